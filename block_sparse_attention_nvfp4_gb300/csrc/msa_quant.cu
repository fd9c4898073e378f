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
// Both roundings equal an exact (real-number) evaluation for every finite input:
//  * scale: the hardware conversion of fl(amax * (1/6)) (relative error below
//    2^-22) is at most one code away from the exact rounding; it is corrected by
//    comparing amax with 6 x the midpoints to its neighbours, 6 v +- 3 x the grid
//    spacing (at most 7 significant bits: exact in FP32).
//  * codes: x / scale correctly rounded to FP32 (reciprocal rounded to nearest, one
//    FMA residual and one FMA correction: Markstein's division), then the hardware
//    round-to-nearest-even conversion to E2M1. The double rounding is harmless: with
//    at most 4 significant bits in the scale, the rounded quotient equals an E2M1
//    midpoint (0.25, 0.75, .. 5) only when x / scale equals it exactly, and lies on
//    the same side of every midpoint as the exact quotient.
//
// Layout: one warp per token; lane = 4 consecutive elements of each of the token's 9
// rows (4 K heads, 4 V heads, the index key), 4 lanes = one 16-element group. All 9
// rows' loads are issued before the token's slot is examined. The 32 group scales of
// the 4 K rows (and of the 4 V rows) are rounded once each, lane 8j + g taking row j's
// group g, and handed back to the group's lanes by shuffles.
#include <cstdint>

#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantCtasPerSm = 3;  // 24 warps x 9 rows x 512 B = 110 KB of loads in flight per SM (80 registers)

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
  const uint32_t e = c >> 3, m = c & 7u;
  const float vc = e4m3_value(c);
  // grid spacing at c: 2^(e-10), 2^-9 for the subnormals; the spacing below c is half
  // of it when c is a power of two above the first binade (m = 0, e >= 2). 6 x the
  // midpoints: 6 vc +- 3 x spacing, at most 7 significant bits: exact.
  const float sp = __uint_as_float((e > 0u ? e + 117u : 118u) << 23);
  const float up = c < 126u ? fmaf(6.f, vc, 3.f * sp) : __int_as_float(0x7f800000);
  const float dn = c > 0u ? fmaf(6.f, vc, (m == 0u && e >= 2u) ? -1.5f * sp : -3.f * sp) : -1.f;
  if (amax > up || (amax == up && (c & 1u))) ++c;
  else if (amax < dn || (amax == dn && (c & 1u))) --c;
  return c;
}

// x / sv correctly rounded, given inv = 1 / sv rounded to nearest; the sign is put back
// for x = -0.0, whose correction step would give +0.0 (-0 + +0 = +0).
__device__ __forceinline__ float div_rn(float x, float sv, float inv) {
  const float q = x * inv;
  return copysignf(fmaf(fmaf(-q, sv, x), inv, q), x);
}

// Two E2M1 codes (sign in bit 3) of x0 / sv (low nibble) and x1 / sv (high nibble).
__device__ __forceinline__ uint32_t e2m1x2(float x0, float x1, float sv, float inv) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r)
      : "f"(div_rn(x1, sv, inv)), "f"(div_rn(x0, sv, inv)));
  return r & 0xFFu;
}

// Largest magnitude of this lane's 16-element group (4 lanes, 4 elements each).
__device__ __forceinline__ float group_amax(const float4& x) {
  float a = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
  return fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
}

// Codes of this lane's 4 elements given its group's scale value and reciprocal, and the
// stores: 2 code bytes per lane, the scale byte by lane 4g.
__device__ __forceinline__ void codes_store(const float4& x, uint32_t sc, float sv, float inv, uint8_t* codes,
                                            uint8_t* scales, int lane) {
  uint32_t c = e2m1x2(x.x, x.y, sv, inv) | (e2m1x2(x.z, x.w, sv, inv) << 8);
  if (sv == 0.f) c = 0u;  // a zero scale gives zero codes
  reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(c);
  if ((lane & 3) == 0) scales[lane >> 2] = static_cast<uint8_t>(sc);
}

// Quantise one 128-element row (this lane's 4 elements) and store it.
__device__ __forceinline__ void quantize_store(const float4& x, uint8_t* codes, uint8_t* scales, int lane) {
  const uint32_t sc = scale_code(group_amax(x));
  const float sv = e4m3_value(sc);
  codes_store(x, sc, sv, __frcp_rn(sv), codes, scales, lane);
}

// Four rows at once: their 32 group scales are rounded once each, lane 8j + g taking
// row j's group g, then handed back to the 4 lanes of each group (the rounding and the
// reciprocal are most of a row's work when every lane repeats them).
__device__ __forceinline__ void quantize_store4(const float4 (&x)[4], uint8_t* const (&codes)[4],
                                                uint8_t* const (&scales)[4], int lane) {
  float am[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) am[j] = group_amax(x[j]);
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float t = __shfl_sync(0xFFFFFFFFu, am[j], 4 * (lane & 7));
    if ((lane >> 3) == j) a = t;
  }
  const uint32_t sc = scale_code(a);
  const float sv = e4m3_value(sc);
  const float inv = __frcp_rn(sv);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int src = 8 * j + (lane >> 2);
    codes_store(x[j], __shfl_sync(0xFFFFFFFFu, sc, src), __shfl_sync(0xFFFFFFFFu, sv, src),
                __shfl_sync(0xFFFFFFFFu, inv, src), codes[j], scales[j], lane);
  }
}

__global__ void __launch_bounds__(kQuantThreads, kQuantCtasPerSm) kv_insert_kernel(const KvInsertParams p) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kQuantThreads / 32);
  for (long long t = static_cast<long long>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
       t < p.num_tokens; t += nwarps) {
    const long long sl = p.slot_mapping[t];
    float4 xk[kGroups], xv[kGroups], xi;
    if (p.k != nullptr)
#pragma unroll
      for (int h = 0; h < kGroups; ++h) xk[h] = __ldcs(reinterpret_cast<const float4*>(p.k + (t * kGroups + h) * kDim) + lane);
    if (p.v != nullptr)
#pragma unroll
      for (int h = 0; h < kGroups; ++h) xv[h] = __ldcs(reinterpret_cast<const float4*>(p.v + (t * kGroups + h) * kDim) + lane);
    if (p.ki != nullptr) xi = __ldcs(reinterpret_cast<const float4*>(p.ki + t * kDim) + lane);
    if (sl < 0) continue;
    const long long page = sl >> 7, slot = sl & 127;
    if (page >= p.num_pages) {
      if (lane == 0) set_flag(p.flags, kFlagBadSlot);
      continue;
    }
    const long long kv_row = page * kGroups * kBlock + slot;  // + h * kBlock for KV head h
    static_assert(kGroups == 4, "the 4 KV heads are quantised together");
    if (p.k != nullptr) {
      uint8_t* const c[4] = {p.k_data + kv_row * 64, p.k_data + (kv_row + kBlock) * 64,
                             p.k_data + (kv_row + 2 * kBlock) * 64, p.k_data + (kv_row + 3 * kBlock) * 64};
      uint8_t* const sc[4] = {p.k_scale + kv_row * 8, p.k_scale + (kv_row + kBlock) * 8,
                              p.k_scale + (kv_row + 2 * kBlock) * 8, p.k_scale + (kv_row + 3 * kBlock) * 8};
      quantize_store4(xk, c, sc, lane);
    }
    if (p.v != nullptr) {
      uint8_t* const c[4] = {p.v_data + kv_row * 64, p.v_data + (kv_row + kBlock) * 64,
                             p.v_data + (kv_row + 2 * kBlock) * 64, p.v_data + (kv_row + 3 * kBlock) * 64};
      uint8_t* const sc[4] = {p.v_scale + kv_row * 8, p.v_scale + (kv_row + kBlock) * 8,
                              p.v_scale + (kv_row + 2 * kBlock) * 8, p.v_scale + (kv_row + 3 * kBlock) * 8};
      quantize_store4(xv, c, sc, lane);
    }
    if (p.ki != nullptr) {
      const long long ki_row = page * kBlock + slot;
      quantize_store(xi, p.ki_data + ki_row * 64, p.ki_scale + ki_row * 8, lane);
    }
  }
}

}  // namespace

cudaError_t launch_kv_insert(const KvInsertParams& prm, int sm_count, cudaStream_t st) {
  const long long blocks_needed = (prm.num_tokens + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  const long long cap = static_cast<long long>(sm_count) * kQuantCtasPerSm;  // one full wave
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  if (grid <= 0) return cudaSuccess;
  kv_insert_kernel<<<grid, kQuantThreads, 0, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace msa
