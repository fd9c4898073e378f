// Device-side building blocks shared by the libmsa kernels: constants, the
// workspace layout, bounded mbarrier waits, TMA / bulk-copy issue, tcgen05
// (TMEM) wrappers, the NVFP4 -> E4M3 dequantisers and the warp top-k.
//
// Sources for the method (cited by tag):
//   [vLLM-zh] vLLM day-0 blog post on MiniMax-M3.1-Flash (Chinese rewrite,
//             agentlenshq.com): "How MiniMax sparse attention works", "Blackwell
//             MSA kernels / dequantising NVFP4 to FP8 with QMUL4", "AMD NVFP4
//             MSA kernel via table lookup".
//   [MSA-fig] "MiniMax goes sparse: reading the M3 attention mechanism from one
//             diagram" (atlascloud.ai), section 1.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

constexpr int kGroups = 4;        // KV heads = GQA groups
constexpr int kHeads = 32;        // query heads
constexpr int kQPerKV = 8;
constexpr int kDim = 128;
constexpr int kBlock = 128;       // tokens per page / KV block
constexpr int kTopK = 16;
constexpr int kMaxRows = 8;       // query rows per request (speculative decode)
constexpr int kMaxReqs = 4096;      // per-request tables live in shared memory

// device error flags (match MSA_FLAG_* in msa.h)
constexpr uint32_t kFlagBadPage = 0x1u;
constexpr uint32_t kFlagBadLength = 0x2u;
constexpr uint32_t kFlagTimeout = 0x4u;
constexpr uint32_t kFlagBadIds = 0x8u;
constexpr uint32_t kFlagBadSlot = 0x10u;

// bounded waits give up after this long (ns of %globaltimer)
constexpr long long kWaitLimitNs = 1000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_flag(uint32_t* flags, uint32_t f) { atomicOr(flags, f); }

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Three-input maximum (one instruction; NaN inputs are ignored as by max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar), "r"(tx)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, for at most kWaitLimitNs.
// On timeout sets the timeout flag and returns false.
static __device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* flags) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = global_ns();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      set_flag(flags, kFlagTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u1(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// Bring [src, src + bytes) into L2 without waiting (bytes a multiple of 16, src 16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits for all of them (release /
// acquire: shared-memory writes before the barrier are visible to the cluster after it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_cluster_u64(uint32_t caddr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(caddr) : "memory");
  return v;
}
__device__ __forceinline__ float ld_cluster_f1(uint32_t caddr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
  return v;
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// Zeros into 16 consecutive TMEM columns of the warp's lanes.
__device__ __forceinline__ void tmem_zero16(uint32_t taddr) {
  const uint32_t z = 0u;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, "
      "%1};" ::"r"(taddr),
      "r"(z)
      : "memory");
}
// tmem_ld32 that also reduces: returns the maximum of this lane's 32 loaded FP32
// columns (NaN ignored, as max.f32 does), computed by the tensor-memory load path
// instead of the ALU. The loaded values themselves are not needed by the callers.
__device__ __forceinline__ float tmem_ld32_max(uint32_t taddr) {
  uint32_t v[32];
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=f"(m)
      : "r"(taddr)
      : "memory");
  return m;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}
// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle. Each K row
// holds 128 bytes of the MN dimension (one swizzle atom); further atoms along MN
// are `mn_atom_bytes` apart (leading byte offset), 8-row K groups 1024 bytes
// apart (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t mn_atom_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((mn_atom_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
// Instruction descriptor, kind::f8f6f4: E4M3 x E4M3 -> F32, K-major A; B K-major
// (b_mn = false: B stored as N rows of K) or MN-major (b_mn = true: K rows of N).
__device__ __forceinline__ uint32_t idesc_e4m3_f32(int M, int N, bool negate_b, bool b_mn = false) {
  return (1u << 4) | (negate_b ? (1u << 14) : 0u) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// D[tmem] (+)= A[tmem] x B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f8_tmemA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p; }" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Weight-stationary form (tcgen05.mma.ws), both operands in shared memory. With
// M = 32 and N = 128 (measured on GB300), D row r is in TMEM lane 32q + r of every
// quadrant q, which holds D columns 32q .. 32q + 31 in 32 TMEM columns from d_tmem.
__device__ __forceinline__ void mma_f8_ws(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.ws.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Weight-stationary form with F16 operands (K = 16 per instruction), both in shared memory.
__device__ __forceinline__ void mma_f16_ws(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.ws.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor, kind::f16: F16 x F16 -> F32, K-major A, B K- or MN-major.
__device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N, bool b_mn) {
  return (1u << 4) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// D[tmem] (+)= A[tmem] x B[smem], F16 operands (K = 16 per instruction).
__device__ __forceinline__ void mma_f16_tmemA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- NVFP4 -> E4M3
// [vLLM-zh, Blackwell kernels] the cache is NVFP4 while queries are FP8, so the
// kernels turn NVFP4 into FP8 before an FP8 MMA. The FP8 value of an element is
// its E2M1 value times its E4M3 group scale, rounded to E4M3. With 256 possible
// scales and 8 E2M1 magnitudes that is a table ([vLLM-zh, AMD NVFP4 MSA kernel
// via table lookup]: 256 scales x 8 magnitudes, pre-rounded to FP8). Here each
// CTA builds it in shared memory with the hardware conversions and byte-permute
// instructions do four lookups at a time.

__device__ __forceinline__ uint32_t cvt_e2m1x2_scaled(uint32_t byte_pair, uint32_t scale_h2) {
  uint32_t h;
  uint16_t e;
  asm("{ .reg .b8 b; cvt.u8.u32 b, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(h) : "r"(byte_pair));
  asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(scale_h2));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e) : "r"(h));
  return e;
}
__device__ __forceinline__ uint32_t e4m3_to_h2_bcast(uint32_t sbyte) {
  uint32_t h;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "r"(sbyte));
  return (h & 0xFFFFu) | (h << 16);
}
// E4M3 images of the magnitudes of E2M1 codes 0..7 times the scale magnitude
// (E4M3 byte s, sign ignored): .x = codes 0..3, .y = codes 4..7, byte k = code k
// (the e2m1x2 conversions take code pairs).
__device__ __forceinline__ uint2 lut_magnitudes(uint32_t s) {
  const uint32_t sc = e4m3_to_h2_bcast(s & 0x7Fu);
  return make_uint2(cvt_e2m1x2_scaled(0x10, sc) | (cvt_e2m1x2_scaled(0x32, sc) << 16),
                    cvt_e2m1x2_scaled(0x54, sc) | (cvt_e2m1x2_scaled(0x76, sc) << 16));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Signed form: 8 elements of code word w (element k in nibble k) -> two words of
// E4M3 bytes, r0 = elements 0..3, r1 = elements 4..7. Magnitudes come from the
// scale's entry (selector bit 3 cleared); the sign of nibble k lands on bit 7 of
// output byte k.
__device__ __forceinline__ void dq8_signed(uint32_t w, uint32_t L0, uint32_t L1, uint32_t& r0, uint32_t& r1) {
  const uint32_t sel = w & 0x77777777u;
  const uint32_t m0 = prmt(L0, L1, sel);
  const uint32_t m1 = prmt(L0, L1, sel >> 16);
  const uint32_t u = w << 4;
  const uint32_t s0 = prmt(w, u, 0x1504);  // byte k's msb = sign of nibble k, k = 0..3
  const uint32_t s1 = prmt(w, u, 0x3726);  // nibbles 4..7
  r0 = m0 ^ (s0 & 0x80808080u);
  r1 = m1 ^ (s1 & 0x80808080u);
}


// ---------------------------------------------------------------- top-k
// [vLLM-zh §How; MSA-fig §1 TopK] One warp selects the blocks of one group:
// the most recent block (nb-1) plus the 15 best of blocks 0..nb-2 by score,
// ties to the lower id; every block when nb <= 16. ids_out gets 16 ascending
// ids, -1 padded. S[c] is block c's score (16-byte aligned rows; plain loads, or
// with kL2 loads that bypass L1 for scores an earlier kernel wrote).
//
// Ranking key: the score's order-preserving integer image in the high word and
// the complemented block id in the low word, so larger key = higher score, then
// lower id; NaN ranks below everything. -0.0 and +0.0 are equal scores (they tie,
// and the lower id wins), so both map to the image of +0.0.
__device__ __forceinline__ uint64_t topk_key(float v, int id) {
  const uint32_t u = v == 0.f ? 0u : __float_as_uint(v);
  uint32_t hi;
  if (v != v) hi = 0u;
  else hi = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(hi) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ int topk_id(uint64_t key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Warp-wide descending bitonic sort of one u64 per lane.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = shfl_xor_u64(v, j);
      const bool up = (lane & k) == 0;          // this k-block sorts descending
      const bool lower = (lane & j) == 0;       // this lane keeps the larger when descending
      const bool keep_max = (up == lower);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// Descending order of a bitonic sequence held one value per lane (half-cleaners only).
__device__ __forceinline__ uint64_t warp_bitonic_merge_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = shfl_xor_u64(v, j);
    const bool lower = (lane & j) == 0;
    v = lower ? (o > v ? o : v) : (o < v ? o : v);
  }
  return v;
}

// The 32 largest of two descending lists (one value per lane), descending: the larger of
// a[i] and b[31 - i] over all i are those 32 values, and they form a bitonic sequence.
__device__ __forceinline__ uint64_t top32_union(uint64_t a, uint64_t b) {
  const int lane = threadIdx.x & 31;
  const uint64_t r = shfl_u64(b, 31 - lane);
  return warp_bitonic_merge_desc(a > r ? a : r);
}

// Keys of candidates c0 .. c1-1 of S (block scores an earlier kernel or another CTA wrote:
// loads bypass L1), id field = candidate index; batch `base` gives lane l the candidates
// c0 + base + 32u + l, u < 8. All 8 loads are issued before the keys are formed.
__device__ __forceinline__ void load_keys8(const float* S, int c0, int c1, int base, uint64_t (&k)[8]) {
  const int lane = threadIdx.x & 31;
  float v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = c0 + base + 32 * u + lane;
    v[u] = c < c1 ? __ldcg(S + c) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = c0 + base + 32 * u + lane;
    k[u] = c < c1 ? topk_key(v[u], c) : 0ull;
  }
}

// Gather the keys >= T of one batch into surv (up to 64), counting all of them.
__device__ __forceinline__ void keep_survivors(const uint64_t (&k)[8], uint64_t T, uint64_t* surv, int& count) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const bool keep = k[u] != 0ull && k[u] >= T;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
    const int pos = count + __popc(bal & ((1u << lane) - 1u));
    if (keep && pos < 64) surv[pos] = k[u];
    count += __popc(bal);
  }
}

// [vLLM-zh §How; MSA-fig §1 TopK] The 15 largest keys of candidates c0 .. c1-1 by one
// warp, descending: lane i < 15 returns the i-th (0 past the end). The 15th largest lane
// maximum T is at most the 15th largest key (the 15 largest lane maxima are 15 distinct
// candidates), so the keys >= T hold the answer; they are gathered (up to 64; scratch
// surv) and sorted. If more than 64 pass (ties), the candidates >= T are merged 32 at a
// time into a running top 32 instead. Ranges of at most 256 candidates are read once,
// into registers; longer ones are streamed twice.
static __device__ __noinline__ uint64_t warp_best15(const float* S, int c0, int c1, uint64_t* surv) {
  constexpr int L = kTopK - 1;
  const int lane = threadIdx.x & 31;
  const int n = c1 - c0;
  uint64_t lmax = 0ull;
  uint64_t kr[8];
  if (n <= 256) {
    load_keys8(S, c0, c1, 0, kr);
#pragma unroll
    for (int u = 0; u < 8; ++u) lmax = kr[u] > lmax ? kr[u] : lmax;
  } else {
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      load_keys8(S, c0, c1, base, k);
#pragma unroll
      for (int u = 0; u < 8; ++u) lmax = k[u] > lmax ? k[u] : lmax;
    }
  }
  const uint64_t T = shfl_u64(warp_sort_desc(lmax), L - 1);
  int count = 0;
  if (n <= 256) {
    keep_survivors(kr, T, surv, count);
  } else {
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      load_keys8(S, c0, c1, base, k);
      keep_survivors(k, T, surv, count);
    }
  }
  __syncwarp();
  uint64_t top;
  if (count <= 32) {
    top = warp_sort_desc(lane < count ? surv[lane] : 0ull);
  } else if (count <= 64) {
    const uint64_t a = warp_sort_desc(surv[lane]);
    const uint64_t b = warp_sort_desc(lane + 32 < count ? surv[lane + 32] : 0ull);
    top = top32_union(a, b);
  } else {
    top = 0ull;
    for (int base = 0; base < n; base += 256) {
      uint64_t k[8];
      if (n <= 256) {
#pragma unroll
        for (int u = 0; u < 8; ++u) k[u] = kr[u];
      } else {
        load_keys8(S, c0, c1, base, k);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t kk = k[u] >= T ? k[u] : 0ull;
        if (__any_sync(0xFFFFFFFFu, kk != 0ull)) top = top32_union(top, warp_sort_desc(kk));
      }
    }
  }
  __syncwarp();
  return lane < L ? top : 0ull;
}

// The 15 best keys of candidates lo .. hi-1 of S by four warps q = 0..3 (128 threads
// meeting at named barrier bar_id): warp q takes a quarter with warp_best15 and warp 0
// merges the four lists (each the exact best 15 of its quarter, so their union holds the
// best 15 of the range). Returns the i-th best key on lane i < 15 of warp 0 (0 past the
// end and on the other warps). Scratch: lists [4][16], surv [4][64].
__device__ __forceinline__ uint64_t quad_best15(const float* S, int lo, int hi, int q, int bar_id, uint64_t* lists,
                                                uint64_t* surv) {
  const int lane = threadIdx.x & 31;
  const int n = hi - lo;
  const int a = lo + q * n / 4, b = lo + (q + 1) * n / 4;
  const uint64_t k = warp_best15(S, a, b, surv + 64 * q);
  if (lane < kTopK) lists[kTopK * q + lane] = k;
  named_bar_sync(bar_id, 128);
  if (q != 0) return 0ull;
  uint64_t top = lane < kTopK ? lists[lane] : 0ull;
#pragma unroll
  for (int w = 1; w < 4; ++w) top = top32_union(top, lane < kTopK ? lists[kTopK * w + lane] : 0ull);
  return lane < kTopK - 1 ? top : 0ull;
}

// The selection of one group from its 15 best candidate keys (one per lane i < 15 of a
// warp, nonzero) and the recent block nb - 1: the 16 ids ascending into ids_out.
__device__ __forceinline__ void write_selection(uint64_t best, int nb, int32_t* ids_out) {
  const int lane = threadIdx.x & 31;
  const int my_id = lane < kTopK - 1 ? topk_id(best) : nb - 1;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    const int other = __shfl_sync(0xFFFFFFFFu, my_id, j);
    rank += other < my_id ? 1 : 0;
  }
  if (lane < kTopK) ids_out[rank] = my_id;
}

// Score loads of the top-k: plain loads (scores in shared memory, or written by
// this CTA), or loads that bypass L1 (scores an earlier kernel wrote).
template <bool kL2>
__device__ __forceinline__ float4 topk_ld4(const float* p) {
  return kL2 ? __ldcg(reinterpret_cast<const float4*>(p)) : *reinterpret_cast<const float4*>(p);
}
template <bool kL2>
__device__ __forceinline__ float topk_ld1(const float* p) {
  return kL2 ? __ldcg(p) : *p;
}

// Exact top-(kTopK-1) of nc candidates by insertion into per-lane sorted lists
// and a 15-round warp merge; the fallback when the threshold filter keeps too many.
template <bool kL2>
static __device__ __noinline__ void topk_by_insertion(const float* S, int nc, int32_t* sel) {
  const int lane = threadIdx.x & 31;
  constexpr int L = kTopK - 1;
  uint64_t list[L];
#pragma unroll
  for (int j = 0; j < L; ++j) list[j] = 0ull;
  for (int c = lane; c < nc; c += 32) {
    const uint64_t key = topk_key(topk_ld1<kL2>(S + c), c);
    if (key > list[L - 1]) {
#pragma unroll
      for (int j = L - 1; j > 0; --j) list[j] = (key > list[j - 1]) ? list[j - 1] : ((key > list[j]) ? key : list[j]);
      list[0] = key > list[0] ? key : list[0];
    }
  }
#pragma unroll 1
  for (int k = 0; k < L; ++k) {
    uint64_t best = list[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = shfl_xor_u64(best, off);
      best = o > best ? o : best;
    }
    if (list[0] == best) {  // keys are unique per block id: exactly one lane
#pragma unroll
      for (int j = 0; j < L - 1; ++j) list[j] = list[j + 1];
      list[L - 1] = 0ull;
    }
    if (lane == 0) sel[k] = topk_id(best);
  }
  __syncwarp();
}

// scratch: 64 u64 per warp (shared memory), for the threshold filter's survivors.
// S may be global or shared memory (callers stage large score rows in shared
// memory, where the passes below do not wait on dependent global round trips).
template <bool kL2 = false>
static __device__ __noinline__ void warp_topk(const float* S, int nb, int32_t* ids_out, uint64_t* scratch) {
  const int lane = threadIdx.x & 31;
  if (nb <= kTopK) {
    if (lane < kTopK) ids_out[lane] = lane < nb ? lane : -1;
    return;
  }
  constexpr int L = kTopK - 1;
  const int nc = nb - 1;  // candidates: every block but the recent one
  int32_t* sel = reinterpret_cast<int32_t*>(scratch + 48);  // 15 winners (kept apart from survivors 0..47)
  // 1. each lane's best key; loads issued 8 at a time (4 blocks per 16-byte load)
  constexpr int kBatch = 32 * 4 * 8;
  uint64_t lmax = 0ull;
  for (int base = 0; base < nc; base += kBatch) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = base + (u * 32 + lane) * 4;
      v[u] = c < nc ? topk_ld4<kL2>(S + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = base + (u * 32 + lane) * 4;
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c + q < nc) {
          const uint64_t k = topk_key(e[q], c + q);
          lmax = k > lmax ? k : lmax;
        }
    }
  }
  // 2. the 15th largest lane maximum bounds the answer: the 15 largest lane maxima
  //    are 15 distinct candidates, so the 15th best candidate is at least that large
  const uint64_t T = shfl_u64(warp_sort_desc(lmax), L - 1);
  // 3. survivors: every candidate with key >= T (contains the exact top 15); the scores
  //    are read again 8 loads at a time (one round trip per 1,024 candidates)
  int count = 0;
  for (int base = 0; base < nc; base += kBatch) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = base + (u * 32 + lane) * 4;
      v[u] = c < nc ? topk_ld4<kL2>(S + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = base + (u * 32 + lane) * 4;
      const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t key = topk_key(e[q], c + q);
        const bool keep = c + q < nc && key >= T;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
        const int pos = count + __popc(bal & ((1u << lane) - 1u));
        if (keep && pos < 48) scratch[pos] = key;  // predicated, no divergent branch
        count += __popc(bal);
      }
    }
  }
  __syncwarp();
  if (count > 48) {
    topk_by_insertion<kL2>(S, nc, sel);
  } else if (count <= 32) {
    // 4. the survivors, one per lane, sorted descending: the top 15 are lanes 0..14
    const uint64_t k = warp_sort_desc(lane < count ? scratch[lane] : 0ull);
    if (lane < L) sel[lane] = topk_id(k);
    __syncwarp();
  } else {
    // 4. exact rank among the survivors
    for (int i = lane; i < count; i += 32) {
      const uint64_t k = scratch[i];
      int rank = 0;
      for (int j = 0; j < count; ++j) rank += scratch[j] > k ? 1 : 0;
      if (rank < L) sel[rank] = topk_id(k);
    }
    __syncwarp();
  }
  // 5. the 15 winners plus the recent block, ascending
  int my_id = lane < L ? sel[lane] : nb - 1;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    const int other = __shfl_sync(0xFFFFFFFFu, my_id, j);
    rank += (other < my_id) ? 1 : 0;
  }
  __syncwarp();
  if (lane < kTopK) ids_out[rank] = my_id;
}

}  // namespace msa
