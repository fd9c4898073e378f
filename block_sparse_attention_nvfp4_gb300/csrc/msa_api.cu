// libmsa C ABI: argument validation, work planning, workspace layout and kernel
// launches for the MSA decode path. The entry points and their contracts are
// declared and documented in include/msa.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/msa.h"
#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr size_t kWsAlign = 256;
size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p *= 2;
  return p;
}

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev & 63];
  if (d.device != dev) {
    int sms = 0, maj = 0, mi = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
    d.sm_count = sms;
    d.major = maj;
    d.minor = mi;
    d.device = dev;
  }
  *out = d;
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

}  // namespace

// 2-D view of an NVFP4 code plane [rows][64 bytes], boxes of 128 rows, 64-byte swizzle.
msa_status encode_code_map(CUtensorMap* map, const uint8_t* base, long long rows) {
  if (get_encode_fn() != cudaSuccess) return MSA_ERR_CUDA;
  cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlock)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_ERR_CUDA;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Host-side checks of everything the host can see. Device-visible values
// (lengths, page ids) are checked by the kernels.
msa_status validate(const msa_decode_args* a, bool need_kv, bool need_idx) {
  if (a == nullptr) return MSA_ERR_INVALID_ARG;
  if (a->num_kv_heads != kGroups || a->q_per_kv != kQPerKV || a->head_dim != kDim || a->block_size != kBlock ||
      a->top_k != kTopK)
    return MSA_ERR_UNSUPPORTED;
  if (a->num_reqs < 0 || a->num_reqs > kMaxReqs || a->total_rows < 0 || a->max_rows_per_req < 1 ||
      a->max_rows_per_req > kMaxRows || a->num_pages < 1 || a->max_pages_per_req < 1)
    return MSA_ERR_INVALID_ARG;
  if (static_cast<long long>(a->total_rows) > static_cast<long long>(a->num_reqs) * a->max_rows_per_req)
    return MSA_ERR_INVALID_ARG;
  if (static_cast<long long>(a->num_pages) * kGroups * kBlock >= (1LL << 31)) return MSA_ERR_UNSUPPORTED;
  if (!(a->sm_scale > 0.f) || !std::isfinite(a->sm_scale)) return MSA_ERR_INVALID_ARG;
  if (a->num_reqs > 0 && (a->context_lens == nullptr || a->q_indptr == nullptr || a->block_table == nullptr))
    return MSA_ERR_INVALID_ARG;
  const bool rows = a->total_rows > 0;
  if (need_idx && ((rows && a->q_idx == nullptr) || a->ki_data == nullptr || a->ki_scale == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (need_kv && ((rows && a->q == nullptr) || a->k_data == nullptr || a->k_scale == nullptr || a->v_data == nullptr ||
                  a->v_scale == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (need_idx && (!aligned16(a->q_idx) || !aligned16(a->ki_data) || !aligned16(a->ki_scale)))
    return MSA_ERR_INVALID_ARG;
  if (need_kv && (!aligned16(a->q) || !aligned16(a->k_data) || !aligned16(a->k_scale) || !aligned16(a->v_data) ||
                  !aligned16(a->v_scale)))
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

msa_status check_device(int* sm_count) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return MSA_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return MSA_ERR_UNSUPPORTED;
  *sm_count = d.sm_count;
  return MSA_OK;
}

namespace {

struct Ws {
  uint32_t* flags;
  float* block_S;
};

msa_status carve(const msa_decode_args* a, void* ws, size_t ws_bytes, Ws* w) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0) return MSA_ERR_WORKSPACE;
  const WsLayout L = ws_layout(a->num_reqs, a->max_pages_per_req);
  if (ws_bytes < L.total) return MSA_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  w->flags = reinterpret_cast<uint32_t*>(base + L.flags);
  w->block_S = reinterpret_cast<float*>(base + L.block_S);
  return MSA_OK;
}

AttnParams attn_params(const msa_decode_args* a, const Ws& w, const Plan& plan, int32_t* ids, uint16_t* out,
                       float* lse) {
  AttnParams p = {};
  p.num_reqs = a->num_reqs;
  p.num_pages = a->num_pages;
  p.max_pages = a->max_pages_per_req;
  p.total_rows = a->total_rows;
  p.context_lens = a->context_lens;
  p.q_indptr = a->q_indptr;
  p.block_table = a->block_table;
  p.block_ids = ids;
  p.q = a->q;
  p.k_data = a->k_data;
  p.k_scale = a->k_scale;
  p.v_data = a->v_data;
  p.v_scale = a->v_scale;
  p.sm_scale_log2 = a->sm_scale * 1.4426950408889634f;
  p.blocks_per_split = plan.blocks_per_split;
  p.splits = plan.splits;
  p.copies = plan.copies;
  p.max_m = kQPerKV * a->max_rows_per_req;
  p.flags = w.flags;
  p.out = out;
  p.lse = lse;
  return p;
}

}  // namespace

int score_stride(int max_pages) { return (max_pages + 3) / 4 * 4; }

Plan make_plan(int num_reqs, int max_rows_per_req, int sm_count) {
  Plan pl;
  // one attention CTA per SM: the fewest blocks per split that fit the (request, group)
  // x split grid into one wave, but at least 2, so a (request, group)'s splits form a
  // cluster of at most 8 CTAs (the portable cluster size) that merges its partials
  const int pairs = num_reqs * kGroups;
  const int target = sm_count > 0 ? sm_count : 1;
  int bps = pairs > 0 ? pow2_ceil((kTopK * pairs + target - 1) / target) : kTopK;
  if (bps < 2) bps = 2;
  if (bps > kTopK) bps = kTopK;
  pl.blocks_per_split = bps;
  pl.splits = kTopK / bps;
  // 4 copies of the <= 32 query rows down the 128-row tile when every request has at most
  // 4 rows (each thread then takes 32 keys of a block), else 2 copies of <= 64 rows
  pl.copies = max_rows_per_req <= 4 ? 4 : 2;
  return pl;
}

WsLayout ws_layout(int num_reqs, int max_pages) {
  WsLayout L;
  size_t off = 0;
  L.flags = off;
  off = align_up(off + 16);
  L.block_S = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(num_reqs) * kGroups * score_stride(max_pages));
  L.total = off;
  return L;
}

msa_status launch_selection(const msa_decode_args* args, int mode, int32_t* ids, float* scores_out, float* tok,
                            long long stride, uint32_t* flags, float* block_S, int sm_count, cudaStream_t st,
                            bool with_topk, int shard, int nshards, uint64_t* dcp_keys) {
  // the scan's shared memory grows with the request count (its page prefix); the exact-score
  // layout leaves room for about 560 requests within the 227 KB a CTA may opt into
  if (select_smem_bytes(args->num_reqs, mode) > 227 * 1024) return MSA_ERR_UNSUPPORTED;
  if (args->num_reqs == 0) return MSA_OK;
  CUtensorMap map;
  msa_status s = encode_code_map(&map, args->ki_data, static_cast<long long>(args->num_pages) * kBlock);
  if (s != MSA_OK) return s;
  SelectParams p = {};
  p.num_reqs = args->num_reqs;
  p.num_pages = args->num_pages;
  p.max_pages = args->max_pages_per_req;
  p.total_rows = args->total_rows;
  p.context_lens = args->context_lens;
  p.q_indptr = args->q_indptr;
  p.block_table = args->block_table;
  p.q_idx = args->q_idx;
  p.ki_scale = args->ki_scale;
  p.block_S = block_S;
  p.s_stride = score_stride(args->max_pages_per_req);
  p.shard = shard;
  p.nshards = nshards;
  p.flags = flags;
  p.block_ids = ids;
  p.block_scores_out = scores_out;
  p.token_scores = tok;
  p.score_stride = stride;
  if (launch_select(map, p, mode, sm_count, st) != cudaSuccess) return MSA_ERR_CUDA;
  if (mode != 1 && with_topk && launch_topk(p, st) != cudaSuccess) return MSA_ERR_CUDA;
  if (dcp_keys != nullptr && launch_dcp_local(p, dcp_keys, st) != cudaSuccess) return MSA_ERR_CUDA;
  return MSA_OK;
}

}  // namespace msa

namespace msa {
namespace {

// One thread waits, through the library's bounded wait, on phase 0 of an mbarrier that
// nothing arrives at: the wait gives up after its limit, sets the timeout flag and returns.
__global__ void selftest_timeout_kernel(uint32_t* flags) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  mbar_fence_init();
  mbar_wait(smem_u32(&bar), 0, flags);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

msa_status msa_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0 || ws_bytes < 256)
    return MSA_ERR_WORKSPACE;
  int sms = 0;
  msa_status s = check_device(&sms);
  if (s != MSA_OK) return s;
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(ws));
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported geometry or device";
    case MSA_ERR_CUDA: return "CUDA runtime error";
    case MSA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MSA_ERR_BAD_TABLE: return "out-of-range page id or length seen on the device";
    case MSA_ERR_TIMEOUT: return "a bounded on-chip wait timed out";
  }
  return "unknown status";
}

msa_status msa_workspace_size(const msa_decode_args* args, size_t* bytes) {
  if (bytes == nullptr) return MSA_ERR_INVALID_ARG;
  msa_status st = validate(args, false, false);
  if (st != MSA_OK) return st;
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return MSA_ERR_CUDA;
  (void)d;
  *bytes = ws_layout(args->num_reqs, args->max_pages_per_req).total;
  return MSA_OK;
}

msa_status msa_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0) return MSA_ERR_WORKSPACE;
  return cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status msa_get_error(void* ws, size_t ws_bytes, void* stream, uint32_t* flags) {
  if (ws == nullptr || ws_bytes < 16 || flags == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
  if (h != 0 && cudaMemsetAsync(ws, 0, sizeof(h), st) != cudaSuccess) return MSA_ERR_CUDA;
  *flags = h;
  if (h & MSA_FLAG_TIMEOUT) return MSA_ERR_TIMEOUT;
  if (h != 0) return MSA_ERR_BAD_TABLE;
  return MSA_OK;
}

static msa_status run_select(const msa_decode_args* args, int mode, int32_t* ids, float* scores_out, float* tok,
                             long long stride, void* ws, size_t ws_bytes, cudaStream_t st) {
  int sms = 0;
  msa_status s = check_device(&sms);
  if (s != MSA_OK) return s;
  if (select_smem_bytes(args->num_reqs, mode) > 227 * 1024) return MSA_ERR_UNSUPPORTED;
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  return launch_selection(args, mode, ids, scores_out, tok, stride, w.flags, w.block_S, sms, st);
}

msa_status msa_index_scores(const msa_decode_args* args, float* scores, int64_t score_stride, void* ws,
                            size_t ws_bytes, void* stream) {
  msa_status s = validate(args, false, true);
  if (s != MSA_OK) return s;
  if (scores == nullptr || score_stride < static_cast<int64_t>(args->max_pages_per_req) * kBlock)
    return MSA_ERR_INVALID_ARG;
  return run_select(args, 1, nullptr, nullptr, scores, score_stride, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

msa_status msa_select_blocks(const msa_decode_args* args, int32_t* block_ids, float* block_scores, void* ws,
                             size_t ws_bytes, void* stream) {
  msa_status s = validate(args, false, true);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr) return MSA_ERR_INVALID_ARG;
  return run_select(args, 0, block_ids, block_scores, nullptr, 0, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

msa_status msa_select_blocks_exact(const msa_decode_args* args, int32_t* block_ids, float* block_scores, void* ws,
                                   size_t ws_bytes, void* stream) {
  msa_status s = validate(args, false, true);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr) return MSA_ERR_INVALID_ARG;
  return run_select(args, 2, block_ids, block_scores, nullptr, 0, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

msa_status msa_dcp_local_topk(const msa_decode_args* args, int32_t rank, int32_t world, uint64_t* cand_keys,
                              void* ws, size_t ws_bytes, void* stream) {
  msa_status s = validate(args, false, true);
  if (s != MSA_OK) return s;
  if (cand_keys == nullptr || (reinterpret_cast<uintptr_t>(cand_keys) & 7u) != 0 || world < 1 ||
      world > MSA_DCP_MAX_WORLD || rank < 0 || rank >= world)
    return MSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((s = check_device(&sms)) != MSA_OK) return s;
  if (select_smem_bytes(args->num_reqs, 0) > 227 * 1024) return MSA_ERR_UNSUPPORTED;
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  return launch_selection(args, 0, nullptr, nullptr, nullptr, 0, w.flags, w.block_S, sms,
                          static_cast<cudaStream_t>(stream), false, rank, world, cand_keys);
}

msa_status msa_dcp_merge_topk(const msa_decode_args* args, int32_t world, int32_t group0, int32_t n_groups,
                              const uint64_t* all_keys, int32_t* block_ids, void* ws, size_t ws_bytes,
                              void* stream) {
  msa_status s = validate(args, false, false);
  if (s != MSA_OK) return s;
  if (all_keys == nullptr || block_ids == nullptr || (reinterpret_cast<uintptr_t>(all_keys) & 7u) != 0 ||
      world < 1 || world > MSA_DCP_MAX_WORLD || group0 < 0 || n_groups < 1 || group0 + n_groups > kGroups)
    return MSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((s = check_device(&sms)) != MSA_OK) return s;
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  if (args->num_reqs == 0) return MSA_OK;
  DcpMergeParams p = {};
  p.num_reqs = args->num_reqs;
  p.max_pages = args->max_pages_per_req;
  p.total_rows = args->total_rows;
  p.context_lens = args->context_lens;
  p.q_indptr = args->q_indptr;
  p.keys = all_keys;
  p.world = world;
  p.group0 = group0;
  p.n_groups = n_groups;
  p.block_ids = block_ids;
  p.flags = w.flags;
  return launch_dcp_merge(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status msa_block_maxpool_topk(const msa_decode_args* args, const float* scores, int64_t score_stride,
                                  int32_t* block_ids, float* block_scores, void* ws, size_t ws_bytes, void* stream) {
  msa_status s = validate(args, false, false);
  if (s != MSA_OK) return s;
  if (scores == nullptr || block_ids == nullptr ||
      score_stride < static_cast<int64_t>(args->max_pages_per_req) * kBlock)
    return MSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((s = check_device(&sms)) != MSA_OK) return s;
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  if (args->num_reqs == 0) return MSA_OK;
  MaxpoolParams p = {};
  p.num_reqs = args->num_reqs;
  p.max_pages = args->max_pages_per_req;
  p.total_rows = args->total_rows;
  p.context_lens = args->context_lens;
  p.q_indptr = args->q_indptr;
  p.scores = scores;
  p.score_stride = score_stride;
  p.block_S = w.block_S;
  p.s_stride = msa::score_stride(args->max_pages_per_req);
  p.block_ids = block_ids;
  p.block_scores_out = block_scores;
  p.flags = w.flags;
  return launch_maxpool_topk(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// fused: the attention kernel selects the ids itself from the block scores the scan left in
// the workspace (and writes them to ids); otherwise it reads the given ids
static msa_status run_attn(const msa_decode_args* args, int32_t* ids, uint16_t* out, float* lse, void* ws,
                           size_t ws_bytes, cudaStream_t st, bool pdl, bool fused, bool small_rows = false) {
  int sms = 0;
  msa_status s = check_device(&sms);
  if (s != MSA_OK) return s;
  const Plan plan = make_plan(args->num_reqs, args->max_rows_per_req, sms);
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  if (args->num_reqs == 0) return MSA_OK;
  // the K and V code planes as [num_pages * 4 * 128 rows][64 bytes] for the tensor copies
  const long long rows = static_cast<long long>(args->num_pages) * kGroups * kBlock;
  CUtensorMap kmap, vmap;
  if ((s = encode_code_map(&kmap, args->k_data, rows)) != MSA_OK) return s;
  if ((s = encode_code_map(&vmap, args->v_data, rows)) != MSA_OK) return s;
  AttnParams p = attn_params(args, w, plan, ids, out, lse);
  if (fused) {
    p.block_S = w.block_S;
    p.s_stride = score_stride(args->max_pages_per_req);
  }
  if (small_rows) return launch_attn_small(kmap, vmap, p, pdl, st) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
  return launch_attn(kmap, vmap, p, pdl, st) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status msa_sparse_attn_decode(const msa_decode_args* args, const int32_t* block_ids, uint16_t* out_bf16,
                                  float* lse, void* ws, size_t ws_bytes, void* stream) {
  msa_status s = validate(args, true, false);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr || out_bf16 == nullptr) return MSA_ERR_INVALID_ARG;
  return run_attn(args, const_cast<int32_t*>(block_ids), out_bf16, lse, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream), false, false);
}

msa_status msa_sparse_attn_decode_small_rows(const msa_decode_args* args, const int32_t* block_ids,
                                             uint16_t* out_bf16, float* lse, void* ws, size_t ws_bytes,
                                             void* stream) {
  msa_status s = validate(args, true, false);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr || out_bf16 == nullptr) return MSA_ERR_INVALID_ARG;
  if (kQPerKV * args->max_rows_per_req > 16) return MSA_ERR_UNSUPPORTED;
  return run_attn(args, const_cast<int32_t*>(block_ids), out_bf16, lse, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream), false, false, true);
}

msa_status msa_decode(const msa_decode_args* args, int32_t* block_ids, uint16_t* out_bf16, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  msa_status s = validate(args, true, true);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr || out_bf16 == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((s = check_device(&sms)) != MSA_OK) return s;
  if (select_smem_bytes(args->num_reqs, 0) > 227 * 1024) return MSA_ERR_UNSUPPORTED;
  Ws w;
  if ((s = carve(args, ws, ws_bytes, &w)) != MSA_OK) return s;
  // the index scan with its block max pool, then the attention, chained by programmatic
  // dependent launch. The top-k runs in a kernel of its own between them (one CTA per
  // request), except (measured on GB300) in two cases where the attention kernel ranks its
  // group's candidates itself, saving a kernel boundary:
  //  * requests may exceed 1,025 blocks and the attention splits each (request, group) over
  //    4 or more CTAs: each CTA of the cluster ranks a share of the candidates and the cluster
  //    merges the shares (one 524,288-token request: 45.5 -> 42-43 us per step);
  //  * every (request, group) is one CTA and no request exceeds 1,025 blocks: the CTA ranks
  //    its group's candidates alone (32 x 65,536 tokens: ~80 -> ~78.5 us per step).
  // Batches with two splits (16 x 131,072) or longer rows in one CTA (64 ragged requests up
  // to 262,144 tokens) are faster with the kernel.
  const Plan plan = make_plan(args->num_reqs, args->max_rows_per_req, sms);
  const bool fused_topk = (args->max_pages_per_req > 1025 && plan.splits >= 4) ||
                          (args->max_pages_per_req <= 1025 && plan.splits == 1);
  if ((s = launch_selection(args, 0, block_ids, nullptr, nullptr, 0, w.flags, w.block_S, sms, st, !fused_topk)) !=
      MSA_OK)
    return s;
  return run_attn(args, block_ids, out_bf16, lse, ws, ws_bytes, st, true, fused_topk);
}

msa_status msa_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t nrows, uint8_t* out_e4m3,
                            int32_t path, void* stream) {
  if (codes == nullptr || scales == nullptr || out_e4m3 == nullptr || nrows < 0 || (path != 0 && path != 1))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 3u) != 0 || (reinterpret_cast<uintptr_t>(out_e4m3) & 3u) != 0)
    return MSA_ERR_INVALID_ARG;
  int sms = 0;
  msa_status s = check_device(&sms);
  if (s != MSA_OK) return s;
  if (nrows == 0) return MSA_OK;
  return launch_dequant_rows(codes, scales, nrows, out_e4m3, path, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}

msa_status msa_kv_insert_nvfp4(const msa_kv_insert_args* a, void* ws, size_t ws_bytes, void* stream) {
  if (a == nullptr || a->num_tokens < 0 || a->num_pages <= 0) return MSA_ERR_INVALID_ARG;
  if (a->num_tokens > 0 && a->slot_mapping == nullptr) return MSA_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if ((a->k != nullptr && (a->k_data == nullptr || a->k_scale == nullptr || misaligned(a->k))) ||
      (a->v != nullptr && (a->v_data == nullptr || a->v_scale == nullptr || misaligned(a->v))) ||
      (a->k_idx != nullptr && (a->ki_data == nullptr || a->ki_scale == nullptr || misaligned(a->k_idx))))
    return MSA_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0 || ws_bytes < kWsAlign)
    return MSA_ERR_WORKSPACE;
  int sms = 0;
  msa_status s = check_device(&sms);
  if (s != MSA_OK) return s;
  if (a->num_tokens == 0 || (a->k == nullptr && a->v == nullptr && a->k_idx == nullptr)) return MSA_OK;
  KvInsertParams p;
  p.num_tokens = a->num_tokens;
  p.num_pages = a->num_pages;
  p.slot_mapping = a->slot_mapping;
  p.k = a->k;
  p.v = a->v;
  p.ki = a->k_idx;
  p.k_data = a->k_data;
  p.k_scale = a->k_scale;
  p.v_data = a->v_data;
  p.v_scale = a->v_scale;
  p.ki_data = a->ki_data;
  p.ki_scale = a->ki_scale;
  p.flags = static_cast<uint32_t*>(ws);
  return launch_kv_insert(p, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
