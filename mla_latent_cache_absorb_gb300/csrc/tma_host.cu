// Host side of the TMA loads: the CUDA driver's tensor-map encoder, looked up once, and the
// encoding of 2D bf16 maps with a small per-thread cache of recent encodings. Kept apart from
// the kernels so that host-only changes leave the kernel sources untouched.
#include "common.cuh"

#include <cudaTypedefs.h>

namespace mla {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once, thread-safely (a function-local static's initialiser runs exactly once)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    if (e != cudaSuccess) (void)cudaGetLastError();   // leave no error of this lookup behind
    return nullptr;
  }();
  return fn;
}

bool make_map_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows, int swizzle_bytes) {
  // The encoding depends only on these arguments, so recent ones are kept per host thread: a
  // decode step encodes up to five maps, mostly the same ones call after call.
  struct Entry {
    const void* base;
    uint64_t inner, rows;
    uint32_t box_inner, box_rows;
    int swizzle;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries];
  thread_local int n_used = 0, next = 0;
  for (int i = 0; i < n_used; ++i) {
    const Entry& en = cache[i];
    if (en.base == base && en.inner == inner && en.rows == rows && en.box_inner == box_inner &&
        en.box_rows == box_rows && en.swizzle == swizzle_bytes) {
      *m = en.map;
      return true;
    }
  }
  if (swizzle_bytes != 128 && swizzle_bytes != 64) return false;
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{base, inner, rows, box_inner, box_rows, swizzle_bytes, *m};
  next = (next + 1) % kEntries;
  if (n_used < kEntries) ++n_used;
  return true;
}

// Rows of C + R bf16 viewed as [rows][C/64 blocks][64]: one box of box_rows rows x box_blocks
// consecutive 64-column blocks lands as box_blocks separate [box_rows][64] tiles, each with the
// 128-byte swizzle (the same image as box_blocks two-dimensional boxes of 64 columns).
bool make_map_row_blocks_bf16(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows,
                              uint32_t n_blocks, uint32_t box_rows, uint32_t box_blocks) {
  struct Entry {
    const void* base;
    uint64_t row_elems, rows;
    uint32_t n_blocks, box_rows, box_blocks;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries];
  thread_local int n_used = 0, next = 0;
  for (int i = 0; i < n_used; ++i) {
    const Entry& en = cache[i];
    if (en.base == base && en.row_elems == row_elems && en.rows == rows && en.n_blocks == n_blocks &&
        en.box_rows == box_rows && en.box_blocks == box_blocks) {
      *m = en.map;
      return true;
    }
  }
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {64, rows, n_blocks};
  cuuint64_t strides[2] = {row_elems * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_blocks};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{base, row_elems, rows, n_blocks, box_rows, box_blocks, *m};
  next = (next + 1) % kEntries;
  if (n_used < kEntries) ++n_used;
  return true;
}

bool tma_encoder_available() { return encode_fn() != nullptr; }

}  // namespace mla
