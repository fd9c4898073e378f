// msa_select_blocks_noalloc: the block selection (index scan with block max
// pool, then top-k) for callers that cannot allocate device memory.
//
// Who needs this: some hosts give a library only the tensors it works on and
// keep the device allocator to themselves (plugin and custom-operator
// interfaces of inference servers, sandboxed extensions), and some decode loops
// must not call cudaMalloc at all, because it can synchronise the device and
// stall every other stream. Such callers cannot provide the workspace that
// msa_select_blocks takes. This entry point runs the same kernels, through the
// same host checks and launch sequence, with their scratch (device error flags,
// block scores) in a fixed buffer compiled into the library instead.
//
// The buffer is kScratchBytes (8 MiB) of device memory that every GPU which
// loads libmsa holds until the process exits. All calls share it, so calls that
// overlap on the GPU (on different streams, or from different host threads)
// race on it and must be serialised by the caller.
#include "../../include/msa.h"
#include "msa_common.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr size_t kFlagsBytes = 256;  // the flags word, padded so the block scores start 256-byte aligned

// The scratch buffer itself. Host code must not use this name as an address:
// it is a host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// Device address of the scratch buffer on the current device. Looked up on every
// call (a lookup, no allocation), so the address stays right if the device's
// context is torn down and made again (cudaDeviceReset), which may move the buffer.
// The first lookup on a device loads the library's device code there if it was not
// loaded yet, which is why the first call on each device should precede any stream
// capture.
cudaError_t scratch_address(uint8_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *out = static_cast<uint8_t*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_select_blocks_noalloc(const msa_decode_args* args, int32_t* block_ids,
                                                float* block_scores, void* stream) {
  msa_status s = validate(args, false, true);
  if (s != MSA_OK) return s;
  if (block_ids == nullptr) return MSA_ERR_INVALID_ARG;
  // scratch layout: error flags (256 B) | block scores [B][4][max_pages rounded up to 4]
  const size_t need = kFlagsBytes + sizeof(float) * static_cast<size_t>(args->num_reqs) * kGroups *
                                        static_cast<size_t>(score_stride(args->max_pages_per_req));
  if (need > kScratchBytes) return MSA_ERR_WORKSPACE;  // the batch needs more than the fixed buffer holds
  int sms = 0;
  if ((s = check_device(&sms)) != MSA_OK) return s;
  uint8_t* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the flags must start at zero (they then report this call's device-side findings);
  // the block maxima are written before they are read
  if (cudaMemsetAsync(base, 0, kFlagsBytes, st) != cudaSuccess) return MSA_ERR_CUDA;
  return launch_selection(args, 0, block_ids, block_scores, nullptr, 0, reinterpret_cast<uint32_t*>(base),
                          reinterpret_cast<float*>(base + kFlagsBytes), sms, st);
}

extern "C" msa_status msa_select_blocks_noalloc_get_error(void* stream, uint32_t* flags) {
  if (flags == nullptr) return MSA_ERR_INVALID_ARG;
  uint8_t* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, base, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
  *flags = h;
  if (h & MSA_FLAG_TIMEOUT) return MSA_ERR_TIMEOUT;
  if (h != 0) return MSA_ERR_BAD_TABLE;
  return MSA_OK;
}
