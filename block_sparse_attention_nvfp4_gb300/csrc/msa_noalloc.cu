// msa_select_blocks_noalloc: the block selection (index scan with block max
// pool, then top-k) for callers that cannot allocate device memory.
//
// Who needs this: some hosts give a library only the tensors it works on and
// keep the device allocator to themselves (plugin and custom-operator
// interfaces of inference servers, sandboxed extensions), and some decode loops
// must not call cudaMalloc at all, because it can synchronise the device and
// stall every other stream. Such callers cannot provide the workspace that
// msa_select_blocks takes. This entry point runs the same kernels with their
// scratch (device error flags, block scores) in a fixed buffer compiled into
// the library instead.
//
// The buffer is kScratchBytes (8 MiB) of device memory that every GPU which
// loads libmsa holds until the process exits. All calls share it, so calls that
// overlap on the GPU (on different streams, or from different host threads)
// race on it and must be serialised by the caller.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/msa.h"
#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;

// The scratch buffer itself. Host code must not use this name as an address:
// it is a host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};  // device address of g_noalloc_scratch, per device

// Device address of the scratch buffer on the current device, looked up once
// per device (the first call on each device does this).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_select_blocks_noalloc(const msa_decode_args* args, int32_t* block_ids,
                                                float* block_scores, void* stream) {
  if (args == nullptr || block_ids == nullptr) return MSA_ERR_INVALID_ARG;
  if (args->num_kv_heads != kGroups || args->q_per_kv != kQPerKV || args->head_dim != kDim ||
      args->block_size != kBlock || args->top_k != kTopK)
    return MSA_ERR_UNSUPPORTED;
  if (args->num_reqs < 0 || args->num_reqs > kMaxReqs || args->total_rows < 0 || args->max_rows_per_req < 1 ||
      args->max_rows_per_req > kMaxRows || args->num_pages < 1 || args->max_pages_per_req < 1 ||
      static_cast<long long>(args->total_rows) > static_cast<long long>(args->num_reqs) * args->max_rows_per_req)
    return MSA_ERR_INVALID_ARG;
  if (static_cast<long long>(args->num_pages) * kGroups * kBlock >= (1LL << 31)) return MSA_ERR_UNSUPPORTED;
  if (args->num_reqs > 0 && (args->context_lens == nullptr || args->q_indptr == nullptr ||
                             args->block_table == nullptr || args->ki_data == nullptr || args->ki_scale == nullptr ||
                             (args->total_rows > 0 && args->q_idx == nullptr)))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(args->q_idx) & 15u) || (reinterpret_cast<uintptr_t>(args->ki_data) & 15u) ||
      (reinterpret_cast<uintptr_t>(args->ki_scale) & 15u))
    return MSA_ERR_INVALID_ARG;

  // scratch layout: error flags (256 B) | block scores [B][4][max_pages rounded up to 4]
  const size_t off_S = 256;
  const size_t need =
      off_S + sizeof(float) * static_cast<size_t>(args->num_reqs) * kGroups * score_stride(args->max_pages_per_req);
  if (need > kScratchBytes) return MSA_ERR_WORKSPACE;  // the batch needs more than the fixed buffer holds

  int dev = 0, maj = 0, mi = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (maj != 10 || mi != 3) return MSA_ERR_UNSUPPORTED;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MSA_ERR_CUDA;
  if (args->num_reqs == 0) return MSA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* s = static_cast<uint8_t*>(base);
  // the flags must start at zero; the block maxima are written before they are read
  if (cudaMemsetAsync(s, 0, off_S, st) != cudaSuccess) return MSA_ERR_CUDA;

  CUtensorMap map;
  {
    // same tensor view of the index-key codes as msa_select_blocks uses
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return MSA_ERR_CUDA;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(args->num_pages) * kBlock};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlock)};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(args->ki_data), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MSA_ERR_CUDA;
  }
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
  p.flags = reinterpret_cast<uint32_t*>(s);
  p.block_S = reinterpret_cast<float*>(s + off_S);
  p.s_stride = score_stride(args->max_pages_per_req);
  p.block_ids = block_ids;
  p.block_scores_out = block_scores;
  if (launch_select(map, p, 0, sms, st) != cudaSuccess) return MSA_ERR_CUDA;
  return launch_topk(p, st) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
