// mla_decode_attn_noalloc: the decode step of mla_decode_attn with its workspace in a fixed
// array of device memory that is part of the library, so the call allocates nothing.
//
// Who needs it: a caller that may not allocate device memory at the moment it decodes. A
// plugin whose host engine owns every byte of device memory and forbids allocation inside
// its execute hook; a server that reserved its whole memory budget at start-up and must not
// grow past it; a latency-bound decode loop that cannot take the device-wide synchronisation
// cudaMalloc/cudaFree imply. Such callers cannot hand mla_decode_attn a workspace sized for
// the batch, so this entry point brings its own.
//
// This is an addition of the library; the descriptions of the method have no counterpart.
#include <cuda_runtime.h>

#include <cstdint>

#include "mla.h"

namespace {

// The whole decode workspace (error word, fused query rows and their residual, split
// partials, merge metadata) lives here. 64 MiB holds, e.g., 128 heads x 64 sequences on a
// 152-SM device; mla_decode_workspace_size says what a given (cfg, B) needs.
__device__ __align__(256) unsigned char g_scratch[MLA_NOALLOC_SCRATCH_BYTES];

// Device address of g_scratch in the current device's context. Looked up on every call, not
// cached: cudaGetSymbolAddress allocates nothing and is cheap once the module is loaded, and
// a cached address would go stale if the context were torn down and recreated (after a
// cudaDeviceReset the module can load at another address).
mla_status scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();   // leave no error behind for the caller's next CUDA call
    return MLA_ERR_CUDA;
  }
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_attn_noalloc(const mla_config* cfg, const void* q, const void* kv_b,
                                              const mla_cache* cache, const int32_t* seq_lens,
                                              const int32_t* positions, float* out, float* lse,
                                              int32_t B, int32_t* device_error, mla_stream_t stream) {
  // size first: a batch the array cannot hold is refused before anything is enqueued
  size_t need = 0;
  mla_status st = mla_decode_workspace_size(cfg, B, &need);
  if (st != MLA_OK) return st;
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  if (device_error != nullptr && (reinterpret_cast<uintptr_t>(device_error) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  void* ws = nullptr;
  st = scratch_address(&ws);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The error word (the first 256 bytes) is the one part of the workspace the kernels read
  // before writing, and it must hold zero when they start: clear it on the stream, every
  // call, so each call reports only its own device errors.
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return MLA_ERR_CUDA;
  st = mla_decode_attn(cfg, q, kv_b, cache, seq_lens, positions, out, lse, B, ws,
                       (size_t)MLA_NOALLOC_SCRATCH_BYTES, stream);
  if (st != MLA_OK) return st;
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
